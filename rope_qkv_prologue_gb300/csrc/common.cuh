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
__device__ __forceinline__ void rope_cos_sin(int32_t pos, uint64_t turns, float* c, float* s) {
  const uint64_t t = static_cast<uint64_t>(static_cast<int64_t>(pos)) * turns;
  const float x = static_cast<float>(static_cast<int64_t>(t)) * 1.0842021724855044e-19f;  // 2^-63
  sincospif(x, s, c);
}

}  // namespace qkvp
