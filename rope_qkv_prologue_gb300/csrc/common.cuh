// Device-side building blocks shared by the prologue kernels (sm_103a).
//
// Data movement: every tensor is moved in 16-byte chunks (8 bf16). A head of
// head_dim = 64 is 8 consecutive chunks, so 8 consecutive lanes of a warp hold
// one head, and the rotate-half partner of element i (element i + D/2) sits in
// lane (lane ^ 4) at the same position of its chunk.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace qkvp {

// -------------------------------------------- programmatic dependent launch ----
//
// Every kernel of the library is launched with programmatic stream
// serialization, so its launch and set-up may overlap the tail of the kernel
// before it in the stream. griddep_wait() blocks until every earlier grid has
// finished and its memory is visible: each kernel calls it before its first
// global-memory access. griddep_launch_dependents() lets the next kernel's
// launch begin (it still waits for this one to finish before touching memory).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::); }

// ---------------------------------------------------------------- bf16 ----

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// --------------------------------------------------------- memory ops ----

// Read-once input stream: cache-streaming load (evict first).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
// Output read soon by the next kernel: plain write-back store.
__device__ __forceinline__ void st_keep(uint4* p, const uint4& v) { *p = v; }
// Output read much later (saved activations): cache-streaming store.
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }

// --------------------------------------------------- paired float math ----
//
// Element-wise math runs on pairs of floats with Blackwell's paired fp32
// instructions (__fmul2_rn / __ffma2_rn: two IEEE float operations, each
// rounded exactly as the scalar operation would be). Every kernel computes a
// chunk through the helpers below, so all code paths (streaming or register,
// contiguous or pool destination) produce the same bits for the same inputs.

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

__device__ __forceinline__ void unpack_pairs(const uint4& v, float2 (&p)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = f2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

__device__ __forceinline__ uint4 pack_pairs(const float2 (&p)[4]) {
  return make_uint4(pack2(p[0].x, p[0].y), pack2(p[1].x, p[1].y), pack2(p[2].x, p[2].y), pack2(p[3].x, p[3].y));
}

__device__ __forceinline__ void load_pairs(const float* p, float2 (&w)[4]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  w[0] = f2(a.x, a.y); w[1] = f2(a.z, a.w); w[2] = f2(b.x, b.y); w[3] = f2(b.z, b.w);
}

// Sum over the CPH lanes of a head of one value per lane, in the head's tree
// order: first each lane with its rotate-half partner (lane ^ CPH/2), then
// xor rounds 1, 2, .., CPH/4. The pair-per-lane kernels hold a chunk and its
// partner in one lane, so they start with a local add and save a round of
// shuffles per sum; the order is the same, so both give the same bits.
template <int CPH>
__device__ __forceinline__ float head_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, CPH / 2);
#pragma unroll
  for (int o = 1; o < CPH / 2; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of squares of this lane's 8 values, then over the CPH lanes of the head.
template <int CPH>
__device__ __forceinline__ float head_sum_sq(const float2 (&x)[4]) {
  float2 a = __fmul2_rn(x[0], x[0]);
  a = __ffma2_rn(x[1], x[1], a);
  a = __ffma2_rn(x[2], x[2], a);
  a = __ffma2_rn(x[3], x[3], a);
  return head_sum<CPH>(a.x + a.y);
}

// x + b on pairs (the qkv bias of the GQAttention variant, added before
// anything else).
__device__ __forceinline__ void add_bias_pairs(float2 (&x)[4], const float2 (&b)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = __fadd2_rn(x[i], b[i]);
}

// Forward of one chunk (8 values of one head, already widened; the head's CPH
// lanes call this together): y = x * r * w with r = (mean(x^2) + eps)^-1/2
// (y = x when NORM is off), then rotate-half: o = y * cos + y_partner * ssin,
// where the partner (element +- D/2) is in lane ^ CPH/2 and ssin = -sin for
// the first half of the head, +sin for the second.
template <int CPH, bool ROPE, bool NORM>
__device__ __forceinline__ void chunk_forward(const float2 (&x)[4], const float2 (&w)[4], float eps, float inv_hd,
                                              const float2 (&c)[4], const float2 (&ssin)[4], float2 (&y)[4]) {
  if (NORM) {
    const float r = rsqrtf(fmaf(head_sum_sq<CPH>(x), inv_hd, eps));
    const float2 rr = f2(r, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = __fmul2_rn(__fmul2_rn(x[i], rr), w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = x[i];
  }
  if (ROPE) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 yp = f2(__shfl_xor_sync(0xffffffffu, y[i].x, CPH / 2),
                           __shfl_xor_sync(0xffffffffu, y[i].y, CPH / 2));
      y[i] = __ffma2_rn(y[i], c[i], __fmul2_rn(yp, ssin[i]));
    }
  }
}

// Backward of one chunk. d: gradient of the roped output; x: the norm's input.
//   g  = R(theta)^T d = d * cos + d_partner * ssin   (ssin = +sin / -sin for
//        the first / second half of the head: the transpose flips the sign)
//   r  = (mean(x^2) + eps)^-1/2
//   dx = r (w g) - x (r^3 / D) sum(x w g)
// Also returns gx = g * x (the weight gradient is gx * r) and r. Without the
// norm dx = g (x, w, gx and r unused).
template <int CPH, bool ROPE, bool NORM>
__device__ __forceinline__ void chunk_backward(const float2 (&d)[4], const float2 (&x)[4], const float2 (&w)[4],
                                               float eps, float inv_hd, const float2 (&c)[4],
                                               const float2 (&ssin)[4], float2 (&dx)[4], float2 (&gx)[4],
                                               float& r_out) {
  float2 g[4], wg[4];
  if (ROPE) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 dp = f2(__shfl_xor_sync(0xffffffffu, d[i].x, CPH / 2),
                           __shfl_xor_sync(0xffffffffu, d[i].y, CPH / 2));
      g[i] = __ffma2_rn(d[i], c[i], __fmul2_rn(dp, ssin[i]));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) g[i] = d[i];
  }
  if (!NORM) {
#pragma unroll
    for (int i = 0; i < 4; ++i) dx[i] = gx[i] = g[i];
    r_out = 0.f;
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) wg[i] = __fmul2_rn(w[i], g[i]);
  float2 sq = __fmul2_rn(x[0], x[0]), dt = __fmul2_rn(x[0], wg[0]);
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    sq = __ffma2_rn(x[i], x[i], sq);
    dt = __ffma2_rn(x[i], wg[i], dt);
  }
  const float ss = head_sum<CPH>(sq.x + sq.y), dot = head_sum<CPH>(dt.x + dt.y);
  const float r = rsqrtf(fmaf(ss, inv_hd, eps));
  const float kx = r * r * r * dot * inv_hd;
  const float2 rr = f2(r, r), nk = f2(-kx, -kx);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dx[i] = __ffma2_rn(x[i], nk, __fmul2_rn(rr, wg[i]));
    gx[i] = __fmul2_rn(g[i], x[i]);
  }
  r_out = r;
}

// ---------------------------------------------- pair-per-lane variants ----
//
// The same arithmetic with a different lane layout: one lane holds chunk e of
// a head ("lo", values 8e .. 8e+7) and its rotate-half partner chunk e + CPH/2
// ("hi"), so CPH/2 lanes share a head. The head sums are added in exactly the
// tree order of head_sum (lo + hi, then xor rounds 1, 2, .. over the CPH/2
// lanes), and the rotation uses the same operations on the same operands, so
// results are bit-identical to chunk_forward / chunk_backward.

__device__ __forceinline__ float chunk_partial_sq(const float2 (&x)[4]) {
  float2 a = __fmul2_rn(x[0], x[0]);
  a = __ffma2_rn(x[1], x[1], a);
  a = __ffma2_rn(x[2], x[2], a);
  a = __ffma2_rn(x[3], x[3], a);
  return a.x + a.y;
}

// Sum over the head of per-chunk partials p_lo, p_hi held by the CPH/2 lanes.
template <int CPH>
__device__ __forceinline__ float pair_head_sum(float lo, float hi) {
  float v = lo + hi;
#pragma unroll
  for (int o = 1; o < CPH / 2; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Forward of a chunk pair (widened, biased): y = x * r * w (y = x without the
// norm), then o_lo = y_lo cos - y_hi sin, o_hi = y_hi cos + y_lo sin (c, sn:
// cos and sin of the lane's 8 frequencies).
template <int CPH, bool ROPE, bool NORM>
__device__ __forceinline__ void pair_forward(const float2 (&lo)[4], const float2 (&hi)[4], const float2 (&wlo)[4],
                                             const float2 (&whi)[4], float eps, float inv_hd, const float2 (&c)[4],
                                             const float2 (&sn)[4], float2 (&ylo)[4], float2 (&yhi)[4]) {
  if (NORM) {
    const float ss = pair_head_sum<CPH>(chunk_partial_sq(lo), chunk_partial_sq(hi));
    const float r = rsqrtf(fmaf(ss, inv_hd, eps));
    const float2 rr = f2(r, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ylo[i] = __fmul2_rn(__fmul2_rn(lo[i], rr), wlo[i]);
      yhi[i] = __fmul2_rn(__fmul2_rn(hi[i], rr), whi[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ylo[i] = lo[i];
      yhi[i] = hi[i];
    }
  }
  if (ROPE) {
    const float2 neg = f2(-1.f, -1.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 ns = __fmul2_rn(sn[i], neg);
      const float2 a = __ffma2_rn(ylo[i], c[i], __fmul2_rn(yhi[i], ns));
      const float2 b = __ffma2_rn(yhi[i], c[i], __fmul2_rn(ylo[i], sn[i]));
      ylo[i] = a;
      yhi[i] = b;
    }
  }
}

// Backward of a chunk pair (see chunk_backward): g_lo = d_lo cos + d_hi sin,
// g_hi = d_hi cos - d_lo sin, then the RMSNorm backward with the head's r
// (x: the norm's input, widened and biased). Without the norm dx = g.
template <int CPH, bool ROPE, bool NORM>
__device__ __forceinline__ void pair_backward(const float2 (&dlo)[4], const float2 (&dhi)[4], const float2 (&xlo)[4],
                                              const float2 (&xhi)[4], const float2 (&wlo)[4], const float2 (&whi)[4],
                                              float eps, float inv_hd, const float2 (&c)[4], const float2 (&sn)[4],
                                              float2 (&dxlo)[4], float2 (&dxhi)[4], float2 (&gxlo)[4],
                                              float2 (&gxhi)[4], float& r_out) {
  float2 glo[4], ghi[4];
  if (ROPE) {
    const float2 neg = f2(-1.f, -1.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 ns = __fmul2_rn(sn[i], neg);
      glo[i] = __ffma2_rn(dlo[i], c[i], __fmul2_rn(dhi[i], sn[i]));
      ghi[i] = __ffma2_rn(dhi[i], c[i], __fmul2_rn(dlo[i], ns));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      glo[i] = dlo[i];
      ghi[i] = dhi[i];
    }
  }
  if (!NORM) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dxlo[i] = gxlo[i] = glo[i];
      dxhi[i] = gxhi[i] = ghi[i];
    }
    r_out = 0.f;
    return;
  }
  float2 wglo[4], wghi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    wglo[i] = __fmul2_rn(wlo[i], glo[i]);
    wghi[i] = __fmul2_rn(whi[i], ghi[i]);
  }
  float2 sql = __fmul2_rn(xlo[0], xlo[0]), sqh = __fmul2_rn(xhi[0], xhi[0]);
  float2 dtl = __fmul2_rn(xlo[0], wglo[0]), dth = __fmul2_rn(xhi[0], wghi[0]);
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    sql = __ffma2_rn(xlo[i], xlo[i], sql);
    sqh = __ffma2_rn(xhi[i], xhi[i], sqh);
    dtl = __ffma2_rn(xlo[i], wglo[i], dtl);
    dth = __ffma2_rn(xhi[i], wghi[i], dth);
  }
  const float ss = pair_head_sum<CPH>(sql.x + sql.y, sqh.x + sqh.y);
  const float dot = pair_head_sum<CPH>(dtl.x + dtl.y, dth.x + dth.y);
  const float r = rsqrtf(fmaf(ss, inv_hd, eps));
  const float kx = r * r * r * dot * inv_hd;
  const float2 rr = f2(r, r), nk = f2(-kx, -kx);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dxlo[i] = __ffma2_rn(xlo[i], nk, __fmul2_rn(rr, wglo[i]));
    dxhi[i] = __ffma2_rn(xhi[i], nk, __fmul2_rn(rr, wghi[i]));
    gxlo[i] = __fmul2_rn(glo[i], xlo[i]);
    gxhi[i] = __fmul2_rn(ghi[i], xhi[i]);
  }
  r_out = r;
}

// ------------------------------------------------------ MLA latent rows ----
//
// Norm part of an MLA latent row: lane l of a warp holds norm chunks l, l + 32,
// ... (NCL of them, zero beyond norm_chunks). Both latent kernels use these,
// so they agree bit for bit.

template <int NCL>
__device__ __forceinline__ float latent_sum_sq(const uint4 (&xr)[NCL], float2 (&x)[NCL][4]) {
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < NCL; ++m) {
    unpack_pairs(xr[m], x[m]);
    ss += chunk_partial_sq(x[m]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return ss;
}

// r = 1 / sqrt(ss / n + eps) for R = 1, 2 or 4 rows at once; s[j] is this
// lane's partial sum of squares of row j, r[j] comes back in every lane.
// The reduction is latent_sum_sq's xor butterfly (partners 16, 8, 4, 2, 1)
// with rows traded instead of copied: at partner 16 a lane keeps the rows of
// its half (h = lane bit 4) and sends the others, at partner 8 (R = 4) it
// keeps one row of the two (g = lane bit 3). Every addition adds the same two
// values as the butterfly does, so each row's sum and r have the bits
// latent_sum_sq gives, with 2 + 1 + 3 shuffles for four rows instead of 20.
template <int R>
__device__ __forceinline__ void latent_rsqrt_rows(const float (&s)[R], float inv_n, float eps, float (&r)[R]) {
  static_assert(R == 1 || R == 2 || R == 4, "1, 2 or 4 rows");
  const int lane = threadIdx.x & 31;
  const bool h = (lane & 16) != 0, g = (lane & 8) != 0;
  float u;
  if constexpr (R == 4) {
    const float t0 = (h ? s[2] : s[0]) + __shfl_xor_sync(0xffffffffu, h ? s[0] : s[2], 16);
    const float t1 = (h ? s[3] : s[1]) + __shfl_xor_sync(0xffffffffu, h ? s[1] : s[3], 16);
    u = (g ? t1 : t0) + __shfl_xor_sync(0xffffffffu, g ? t0 : t1, 8);  // row 2h + g
  } else if constexpr (R == 2) {
    u = (h ? s[1] : s[0]) + __shfl_xor_sync(0xffffffffu, h ? s[0] : s[1], 16);  // row h
    u += __shfl_xor_sync(0xffffffffu, u, 8);
  } else {
    u = s[0] + __shfl_xor_sync(0xffffffffu, s[0], 16);
    u += __shfl_xor_sync(0xffffffffu, u, 8);
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
  const float rr = rsqrtf(fmaf(u, inv_n, eps));
#pragma unroll
  for (int j = 0; j < R; ++j) r[j] = R == 1 ? rr : __shfl_sync(0xffffffffu, rr, j * (32 / R));
}

__device__ __forceinline__ uint4 latent_norm_chunk(const float2 (&x)[4], float r, const float2 (&w)[4]) {
  const float2 rr = f2(r, r);
  float2 y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = __fmul2_rn(__fmul2_rn(x[i], rr), w[i]);
  return pack_pairs(y);
}

// Rotate-half of one rope chunk pair: lo = values 8e .. 8e+7 of the rope
// part, hi = their partners 8e + 32 .. (c, sn: cos / sin of frequencies
// 8e .. 8e+7).
__device__ __forceinline__ void latent_rope_pair(const uint4& rlo, const uint4& rhi, const float (&c)[8],
                                                 const float (&sn)[8], uint4& olo, uint4& ohi) {
  float xl[8], xh[8], yl[8], yh[8];
  unpack8(rlo, xl);
  unpack8(rhi, xh);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    yl[i] = fmaf(xl[i], c[i], xh[i] * -sn[i]);
    yh[i] = fmaf(xh[i], c[i], xl[i] * sn[i]);
  }
  olo = pack8(yl);
  ohi = pack8(yh);
}

// The same rotation for half a chunk pair: lo = values 8e + 4h .. 8e + 4h + 3
// of the rope part, hi = their partners 32 further on (c, sn: cos / sin of
// those four frequencies).
__device__ __forceinline__ void latent_rope_quad(const uint2& rlo, const uint2& rhi, const float (&c)[4],
                                                 const float (&sn)[4], uint2& olo, uint2& ohi) {
  const float xl[4] = {__uint_as_float(rlo.x << 16), __uint_as_float(rlo.x & 0xffff0000u),
                       __uint_as_float(rlo.y << 16), __uint_as_float(rlo.y & 0xffff0000u)};
  const float xh[4] = {__uint_as_float(rhi.x << 16), __uint_as_float(rhi.x & 0xffff0000u),
                       __uint_as_float(rhi.y << 16), __uint_as_float(rhi.y & 0xffff0000u)};
  float yl[4], yh[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    yl[i] = fmaf(xl[i], c[i], xh[i] * -sn[i]);
    yh[i] = fmaf(xh[i], c[i], xl[i] * sn[i]);
  }
  olo = make_uint2(pack2(yl[0], yl[1]), pack2(yl[2], yl[3]));
  ohi = make_uint2(pack2(yh[0], yh[1]), pack2(yh[2], yh[3]));
}

// ---------------------------------------------------------- division ----

// n / d for n < 2^16 and 2 <= d <= 2^16 with m = floor(2^32 / d) + 1:
// n * m / 2^32 = n / d + n * delta / 2^32 with 0 < delta <= 1, and the error
// term is below 2^-16 <= 1/d, so it never crosses the next integer.
__device__ __forceinline__ uint32_t small_div(uint32_t n, uint32_t m) { return __umulhi(n, m); }

// --------------------------------------------------------------- RoPE ----

// cos and sin of the angle pos * inv_freq, where the angle per unit position
// is held as an unsigned 0.64 fixed-point fraction of a turn
// (turns = frac(inv_freq / 2pi) * 2^64). The product pos * turns modulo 2^64
// is the angle reduced exactly to one turn; read as a signed number it is
// the angle / pi scaled by 2^63, in [-1, 1).
// Both are then multiplied by `scale` (the cos/sin factor of YaRN-style
// scalings; exactly 1 for plain RoPE, which leaves the values unchanged).
__device__ __forceinline__ void rope_cos_sin(int32_t pos, uint64_t turns, float scale, float* c, float* s) {
  const uint64_t t = static_cast<uint64_t>(static_cast<int64_t>(pos)) * turns;
  const float x = static_cast<float>(static_cast<int64_t>(t)) * 1.0842021724855044e-19f;  // 2^-63
  sincospif(x, s, c);
  *c *= scale;
  *s *= scale;
}

}  // namespace qkvp
