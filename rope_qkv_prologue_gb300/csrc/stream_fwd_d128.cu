// Streaming forward kernel instances for head_dim 128.
#include "gqa_stream.cuh"

namespace qkvp {

namespace {
template <bool S, bool R, bool SV, bool P>
const void* ptr() {
  constexpr StreamShape sh = fwd_stream_shape(SV);
  return reinterpret_cast<const void*>(&qkvp_fwd_stream_kernel<128, S, R, SV, P, sh.warps, sh.ctas_per_sm>);
}
template <bool S, bool R>
const void* pick(const FwdVariant& v) {
  if (v.pool) return ptr<S, R, false, true>();
  return v.save_pre ? ptr<S, R, true, false>() : ptr<S, R, false, false>();
}
}  // namespace

const void* fwd_stream_kernel_d128(const FwdVariant& v) {
  if (v.sectioned) return v.rope ? pick<true, true>(v) : pick<true, false>(v);
  return v.rope ? pick<false, true>(v) : pick<false, false>(v);
}

}  // namespace qkvp
